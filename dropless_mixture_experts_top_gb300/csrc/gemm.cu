// gemm.cu -- persistent grouped GEMMs over ragged expert segments on the
// 5th-generation tensor core (tcgen05, sm_103a), one CTA pair per tile.
//
// A grouped GEMM handles every expert's matrix product in one launch, each at
// its real token count, computing only the valid regions; counts stay on the
// device so nothing is copied to the host (NVIDIA MoE article,
// "Optimizacion 1, el GEMM agrupado").  Two shapes of raggedness occur:
//   ragged M  (forward GEMMs, dA, dX): rows = the expert's permuted rows;
//             output tiles of 256 rows start at each expert's first row, rows
//             past the expert's end are computed but never stored.
//   ragged K  (weight gradients): the reduction runs over the expert's rows;
//             each expert gets its own tensor maps whose row extent ends at the
//             expert's last row, so the last 64-row K block is zero-filled past
//             it by the TMA unit itself; an expert with no rows gets an
//             all-zero gradient.
//
// Kernel structure: clusters of two CTAs (a CTA pair on two SMs), persistent,
// static round-robin over 256x256 output tiles.  Each CTA holds 128 rows of A
// and 128 columns of B in a shared-memory ring (3 stages of 128 of K; dA: 5
// stages of 64 of K, its shared memory also holding a G/U ring), so each SM
// reads half the B operand it would need alone; the pair's MMAs (cta_group::2,
// M=256, N=256, K=16, bf16 in, fp32 accumulate) are issued by the first CTA and
// write each CTA's 128 accumulator rows into its own TMEM.
//   warp 0      TMA producer (both CTAs): 128B-swizzled boxes into its ring;
//               both CTAs' copies complete on CTA 0's barrier
//   warp 1      CTA 0: MMA issuer (CTA 1's warp 1 only shares the TMEM allocation)
//   warps 2..    epilogue (both CTAs): tcgen05.ld of its 128 rows from two
//               double-buffered 256-column accumulators, fused SwiGLU /
//               dSwiGLU, bf16 stores; 4 warps (one per TMEM lane quarter), 8
//               (two per quarter, one per column half) for the modes with the
//               heaviest epilogues: gate/up, dA and the router's dx
//   dA only     one more warp streams each tile's G and U into the G/U ring
//   forward GEMMs of an MXFP8 backward: after each tile's epilogue, the
//               epilogue warps quantise part of the weights into the backward's
//               weight codes (8 epilogue warps for the down GEMM too)
// Every wait is bounded; on a timeout the kernel flags the status word,
// drains its own copies and MMAs, frees TMEM and returns.
#include <cuda.h>

#include "common.cuh"
#include "epilogue.cuh"

namespace moe {
namespace {

constexpr int BM = 128;   // rows per CTA (TMEM lanes); a tile is 2*BM rows
constexpr int BN = 256;   // tile columns (TMEM columns per accumulator); BN/2 per CTA
constexpr int BK = 64;    // K per operand box: one 128-byte swizzle row of bf16
constexpr int kABox = BM * BK * 2;            // 16 KB: this CTA's rows of A for 64 of K
constexpr int kBBox = (BN / 2) * BK * 2;      // 16 KB: this CTA's columns of B for 64 of K
// A pipeline stage holds HALVES consecutive 64-wide K blocks of both operands
// ([A k0 | A k1 | B k0 | B k1]): 128 of K, so eight MMAs per barrier round
// trip; dA keeps 64 (its shared memory also holds the G/U ring).
__host__ __device__ constexpr int halves_of(int mode) { return mode == kBwdDA ? 1 : 2; }
__host__ __device__ constexpr int stage_bytes(int mode) { return halves_of(mode) * (kABox + kBBox); }
constexpr int kBox = 64 * 64 * 2;             // one 64x64 bf16 box (MN-major pieces)
constexpr int kMapsPerExpert = 3;             // ragged K: A, B0, B1
// Warps: producer, MMA issuer, then 4 epilogue warps (one per TMEM lane
// quarter).  The epilogue-heavy modes run 8 (two per quarter, one per column
// half): gate/up writes four outputs per element, dA's dSwiGLU reads G and U
// and writes dG and dU, and the router's dx reads and rewrites dx after a
// K = E reduction too short to hide it -- dA also has a warp that streams each
// tile's G and U into a shared-memory ring ahead of its epilogue, and an
// operand ring of 5 stages to make room.  The other modes run slower with 8
// epilogue warps.
__host__ __device__ constexpr int stages_of(int mode) { return mode == kBwdDA ? 5 : 3; }
__host__ __device__ constexpr int epi_warps(int mode, bool wq = false) {
  return (mode == kBwdDA || mode == kFwdGateUp || mode == kRouterDX || (mode == kFwdDown && wq)) ? 8 : 4;
}
__host__ __device__ constexpr int gu_warps(int mode) { return mode == kBwdDA ? 1 : 0; }
__host__ __device__ constexpr int threads_of(int mode, bool wq = false) {
  return 64 + 32 * (epi_warps(mode, wq) + gu_warps(mode));
}
constexpr uint32_t kTmemCols = 2 * BN;
// Shared memory (from a 1024-aligned base): operand stages | barriers (512) |
// three [E+1] tables | epilogue staging tiles | dA: the G/U ring (1024-aligned).
__host__ __device__ constexpr int epi_off(int mode) {
  return (stages_of(mode) * stage_bytes(mode) + 512 + 3 * (kMaxExperts + 1) * 4 + 15) / 16 * 16;
}
__host__ __device__ constexpr int gu_off(int mode, bool wq = false) {
  return (epi_off(mode) + epi_warps(mode, wq) * kEpiTileBytes + 1023) / 1024 * 1024;
}
__host__ __device__ constexpr int smem_bytes(int mode, bool wq = false) {
  return gu_off(mode, wq) + gu_warps(mode) * kGuSlots * kGuChunkBytes + 1024 /*align*/;
}
static_assert(smem_bytes(kBwdDA) <= 227 * 1024 && smem_bytes(kFwdGateUp) <= 227 * 1024 &&
                  smem_bytes(kFwdDown, true) <= 227 * 1024,
              "shared memory budget");

struct Params {
  int M_rows, H, I, E;
  const int32_t *offsets;
  const uint16_t *G, *U;  // dSwiGLU epilogue inputs
  const float *w_row;     // router weight of each permuted row
  float *g_part;          // dA: partial router-weight gradients [M][g_np] (or null)
  int g_np;               // dA: partials per row (2 per 256-column tile)
  uint16_t *o0, *o1, *o2, *o3;
  uint8_t *aw_t, *aw_t_sf;  // gate/up for an MXFP8 backward: w * A along tokens [I, Mpad] (or null)
  int Mpad;
  // forward GEMMs for an MXFP8 backward: the bf16 weights ([E*H, I] gate (0) and
  // up (1), or [E*I, H] down (0)) and their codes along the last axis with scale atoms
  const uint16_t *wsrc[2];
  uint8_t *wq[2], *wq_sf[2];
  float *of;   // router projection: fp32 output
  int n_out;   // router projection: output columns (E)
  int32_t *status;
  const CUtensorMap *expert_maps;  // ragged K: [E][kMapsPerExpert] maps ending at each expert's end
  int kdim;     // ragged M: the fixed reduction length
  int n_tiles;  // column tiles per row tile
  int m_tiles;  // ragged K: row tiles per expert
};

template <int MODE>
struct Traits {
  static constexpr bool kRaggedK = (MODE == kBwdDWDown || MODE == kBwdDWGateUp || MODE == kRouterDW);
  static constexpr int kAMN = kRaggedK ? 1 : 0;  // A operand MN-major in smem
  static constexpr int kBMN =
      (MODE == kFwdGateUp || MODE == kFwdDown || MODE == kRouterFwd || kRaggedK) ? 1 : 0;
  // column tile = [first source | second source], 128 columns each (gate | up):
  // CTA 0 holds the first source's columns, CTA 1 the second's
  static constexpr bool kPair = (MODE == kFwdGateUp || MODE == kBwdDWGateUp);

  static constexpr uint32_t kIdesc = idesc_bf16(2 * BM, BN, kAMN, kBMN);
};

template <int MODE>
__device__ __forceinline__ Tile decode_tile(int tile, const Params &p, const int *s_tp,
                                            const int *s_off, const int *s_pad) {
  using Tr = Traits<MODE>;
  Tile t;
  if constexpr (!Tr::kRaggedK) {
    const int mt_lin = tile / p.n_tiles, nt = tile % p.n_tiles;
    int lo = 0, hi = p.E - 1;  // largest e with s_tp[e] <= mt_lin
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_tp[mid] <= mt_lin)
        lo = mid;
      else
        hi = mid - 1;
    }
    t.e = lo;
    t.m0 = s_off[lo] + (mt_lin - s_tp[lo]) * (2 * BM);
    t.row_end = s_off[lo + 1];
    t.n0 = nt * (Tr::kPair ? BN / 2 : BN);
    t.nkb = p.kdim / BK;
    // the padded token axis of an MXFP8 backward (each expert from a multiple of 128)
    t.krow0 = s_pad[lo] + (t.m0 - s_off[lo]);
    t.kcount = s_pad[lo] + (s_off[lo + 1] - s_off[lo] + 127) / 128 * 128;
  } else {
    const int per = p.m_tiles * p.n_tiles;
    t.e = s_tp[tile / per];  // experts in decreasing order of rows
    const int rem = tile % per;
    t.m0 = (rem / p.n_tiles) * (2 * BM);
    t.n0 = (rem % p.n_tiles) * (Tr::kPair ? BN / 2 : BN);
    t.krow0 = s_off[t.e];
    t.kcount = s_off[t.e + 1] - s_off[t.e];
    t.nkb = (t.kcount + BK - 1) / BK;
    t.row_end = 0;
  }
  return t;
}

// One box into this CTA's stage, completing on CTA 0's barrier for the stage.
struct StageLoad {
  uint32_t bar_cl;  // CTA 0's full barrier for the stage (shared::cluster address)
  __device__ __forceinline__ void operator()(void *dst, const CUtensorMap *m, int c0, int c1) const {
    tma_load_2d_pair(dst, m, bar_cl, c0, c1);
  }
};

// This CTA's share of one stage: 128 rows of A, 128 columns of B.
// This CTA's rows of A in a ragged M tile: all 128 (one box), or, where the
// expert's rows end inside them, the 32-row boxes that hold its rows (nbox of
// them; the MMA reads the rest of the slot, whose rows are never stored).
template <class Load>
__device__ __forceinline__ void load_a_rows(const Load &ld, uint8_t *sa, const CUtensorMap *full,
                                            const CUtensorMap *part, int k0, int arow, int nbox) {
  if (nbox >= 4) {
    ld(sa, full, k0, arow);
  } else {
    for (int b = 0; b < nbox; ++b) ld(sa + b * 32 * BK * 2, part, k0, arow + 32 * b);
  }
}
__device__ __forceinline__ int a_boxes(const Tile &t, int rank) {
  const int valid = t.row_end - (t.m0 + BM * rank);
  return valid >= BM ? 4 : (valid > 0 ? (valid + 31) / 32 : 0);
}

template <int MODE, class Load>
__device__ __forceinline__ void produce_stage(const Tile &t, int kb, int rank, uint8_t *sa,
                                              uint8_t *sb, const Load &ld, const Params &p,
                                              const CUtensorMap *a0, const CUtensorMap *a1,
                                              const CUtensorMap *b0, const CUtensorMap *b1,
                                              const CUtensorMap *a0s, const CUtensorMap *a1s) {
  const int arow = t.m0 + BM * rank;        // ragged M: this CTA's rows of A
  const int nbox = a_boxes(t, rank);
  const int bcol = t.n0 + (BN / 2) * rank;  // this CTA's columns of B (unpaired modes)
  if constexpr (MODE == kFwdGateUp) {
    load_a_rows(ld, sa, a0, a0s, kb * BK, arow, nbox);
    const CUtensorMap *w = rank == 0 ? b0 : b1;  // gate columns | up columns
    const int wrow = t.e * p.H + kb * BK;
    ld(sb, w, t.n0, wrow);
    ld(sb + kBox, w, t.n0 + 64, wrow);
  } else if constexpr (MODE == kFwdDown || MODE == kRouterFwd) {
    load_a_rows(ld, sa, a0, a0s, kb * BK, arow, nbox);
    const int wrow = t.e * p.I + kb * BK;
    ld(sb, b0, bcol, wrow);
    ld(sb + kBox, b0, bcol + 64, wrow);
  } else if constexpr (MODE == kBwdDA || MODE == kRouterDX) {
    load_a_rows(ld, sa, a0, a0s, kb * BK, arow, nbox);
    ld(sb, b0, kb * BK, t.e * p.I + bcol);
  } else if constexpr (MODE == kBwdDX) {
    const int kbi = p.I / BK;
    if (kb < kbi) {
      load_a_rows(ld, sa, a0, a0s, kb * BK, arow, nbox);
      ld(sb, b0, kb * BK, t.e * p.H + bcol);
    } else {
      load_a_rows(ld, sa, a1, a1s, (kb - kbi) * BK, arow, nbox);
      ld(sb, b1, (kb - kbi) * BK, t.e * p.H + bcol);
    }
  } else if constexpr (MODE == kBwdDWDown || MODE == kRouterDW) {
    const CUtensorMap *em = p.expert_maps + t.e * kMapsPerExpert;  // rows end at the expert's end
    const int r = t.krow0 + kb * BK;
    ld(sa, em + 0, t.m0 + BM * rank, r);
    ld(sa + kBox, em + 0, t.m0 + BM * rank + 64, r);
    ld(sb, em + 1, bcol, r);
    ld(sb + kBox, em + 1, bcol + 64, r);
  } else {  // kBwdDWGateUp
    const CUtensorMap *em = p.expert_maps + t.e * kMapsPerExpert;
    const int r = t.krow0 + kb * BK;
    ld(sa, em + 0, t.m0 + BM * rank, r);
    ld(sa + kBox, em + 0, t.m0 + BM * rank + 64, r);
    const CUtensorMap *g = em + (rank == 0 ? 1 : 2);  // dG columns | dU columns
    ld(sb, g, t.n0, r);
    ld(sb + kBox, g, t.n0 + 64, r);
  }
}

// The backward's weight codes for 32 rows x 128 columns of a bf16 weight
// ([rows, ld] row-major, row0 a multiple of 32, col0 of 128): E4M3 codes and
// UE8M0 scales in blocks of 32 along the rows, the quantiser's rule
// (mxfp8.cuh).  One warp: four rows per step, eight lanes per row, sixteen
// columns per lane, so a block's amax takes one exchange between lane pairs and
// each row leaves as one 128-byte line of codes and one 4-byte word of scales.
// The 32 rows lie in one 128-row scale atom (segments and groups are multiples
// of 64 rows), so the scale words are the atom's base plus the row's offset.
// Each batch of kBatch steps issues its loads together (all eight where the
// kernel's registers allow).
template <int kBatch>
__device__ __forceinline__ void quant_weight_rows(const uint16_t *__restrict__ w, int row0, int col0, int ld,
                                                  uint8_t *__restrict__ codes, uint8_t *__restrict__ sf,
                                                  SfLayout L, int lane) {
  const int sub = lane & 7, r4 = lane >> 3;
  const size_t base = atom_byte(row0, col0 >> 5, ld, L);  // word of the block's first row
  const int w0 = (row0 - (row0 / L.seg) * L.seg) % L.group & 127;  // its row within the atom
  const uint4 *src = reinterpret_cast<const uint4 *>(w + static_cast<size_t>(row0 + r4) * ld + col0 + sub * 16);
  uint8_t *dst = codes + static_cast<size_t>(row0 + r4) * ld + col0 + sub * 16;
  const size_t step = static_cast<size_t>(4) * ld;  // four rows, in elements and in code bytes
#pragma unroll 1
  for (int bt = 0; bt < 8 / kBatch; ++bt) {
    uint4 in[kBatch][2];
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const size_t off = (bt * kBatch + j) * step / 8;
      in[j][0] = __ldg(src + off);
      in[j][1] = __ldg(src + off + 1);
    }
#pragma unroll
    for (int j = 0; j < kBatch; ++j) {
      const int i = bt * kBatch + j;  // step: rows 4i .. 4i+3 of the 32
      const uint32_t u[8] = {in[j][0].x, in[j][0].y, in[j][0].z, in[j][0].w,
                             in[j][1].x, in[j][1].y, in[j][1].z, in[j][1].w};
      float v[16];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        v[2 * q] = bf16_lo(u[q]);
        v[2 * q + 1] = bf16_hi(u[q]);
      }
      float m[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        m[q] = fmaxf(fmaxf(fabsf(v[q]), fabsf(v[q + 4])), fmaxf(fabsf(v[q + 8]), fabsf(v[q + 12])));
      float amax = fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));  // the other half of the block
      const int X = mx_scale_exp(amax);
      const float sc = pow2_neg(X);
      uint4 o;
      o.x = pack_e4m3x4_scaled(v[0], v[1], v[2], v[3], sc);
      o.y = pack_e4m3x4_scaled(v[4], v[5], v[6], v[7], sc);
      o.z = pack_e4m3x4_scaled(v[8], v[9], v[10], v[11], sc);
      o.w = pack_e4m3x4_scaled(v[12], v[13], v[14], v[15], sc);
      *reinterpret_cast<uint4 *>(dst + i * step) = o;
      // the row's four blocks: scale codes of lanes 0, 2, 4, 6 of its eight, one word
      const uint32_t x0 = static_cast<uint32_t>(X + 127);
      const uint32_t x1 = __shfl_down_sync(0xffffffffu, x0, 2);
      const uint32_t x2 = __shfl_down_sync(0xffffffffu, x0, 4);
      const uint32_t x3 = __shfl_down_sync(0xffffffffu, x0, 6);
      if (sub == 0) {
        const int wr = w0 + 4 * i + r4;  // the row within its atom
        *reinterpret_cast<uint32_t *>(sf + base + (wr & 31) * 16 + (wr >> 5) * 4 - (w0 & 31) * 16 - (w0 >> 5) * 4) =
            x0 | (x1 << 8) | (x2 << 16) | (x3 << 24);
      }
    }
  }
}

template <int MODE, bool WQ>
__global__ void __launch_bounds__(threads_of(MODE, WQ), 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA0,
                        const __grid_constant__ CUtensorMap tmA1,
                        const __grid_constant__ CUtensorMap tmB0,
                        const __grid_constant__ CUtensorMap tmB1,
                        const __grid_constant__ CUtensorMap tmA0s,
                        const __grid_constant__ CUtensorMap tmA1s, const Params p) {
  using Tr = Traits<MODE>;
  static_assert(!WQ || MODE == kFwdGateUp || MODE == kFwdDown, "weight codes come from the forward GEMMs");
  constexpr int STAGES = stages_of(MODE), HALVES = halves_of(MODE);
  constexpr int NT = threads_of(MODE, WQ), EW = epi_warps(MODE, WQ);
  constexpr int kStageBytes = stage_bytes(MODE), kABytes = HALVES * kABox;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *stages = smem;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGES * kStageBytes);
  uint64_t *full = bars;                 // [STAGES] CTA 0 only: both CTAs' copies landed
  uint64_t *empty = bars + STAGES;       // [STAGES] pair MMA (and weight quantisers) done with the stage
  uint64_t *tfull = bars + 2 * STAGES;   // [2] accumulator ready (both CTAs)
  uint64_t *tempty = tfull + 2;          // [2] CTA 0 only: both CTAs' epilogues done
  uint64_t *drain = tempty + 2;          // abort path: MMA completion
  uint64_t *gu_full = drain + 1;         // [kGuSlots] dA: a G/U chunk landed (this CTA)
  uint64_t *gu_empty = gu_full + kGuSlots;  // [kGuSlots] dA: its 4 epilogue warps read it
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gu_empty + kGuSlots);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  // [E+1] ragged M: tile prefix over experts; ragged K: experts by decreasing row count
  int *s_tp = reinterpret_cast<int *>(smem + STAGES * kStageBytes + 512);
  int *s_off = s_tp + (kMaxExperts + 1);                                    // [E+1] row offsets
  int *s_pad = s_off + (kMaxExperts + 1);  // [E+1] ragged M: padded offsets (128-aligned segments)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;
  const int rank = static_cast<int>(cluster_ctarank());  // 0: issues the pair's MMAs
  uint8_t *epi_tiles = smem + epi_off(MODE);  // [epilogue warp] 32 x 32 bf16 staging tiles
  uint8_t *gu_ring = smem + gu_off(MODE, WQ); // dA: [kGuSlots] G chunk | U chunk
  const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 2 * EW);  // one arrival per epilogue warp of both CTAs
    }
    mbar_init(drain, 1);
    for (int s = 0; s < kGuSlots; ++s) {
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
  if (warp == 1) tmem_alloc_pair(tmem_slot, kTmemCols);
  griddep_wait();  // the set-up above overlaps the previous kernel's end; its outputs are read below
  // no offsets: one segment of all M_rows rows (the router projection's logits and dx)
  for (int e = threadIdx.x; e <= E; e += NT)
    s_off[e] = p.offsets ? __ldg(p.offsets + e) : (e == 0 ? 0 : p.M_rows);
  __syncthreads();
  bool skewed = false;
  if (Tr::kRaggedK) {
    // Skewed routing (an expert with more than twice the mean rows): longest
    // reductions first, and the tiles go out in a snake over the CTA pairs
    // (round r to pairs 0, 1, ... when r is even, to pairs ..., 1, 0 when odd),
    // which balances decreasing work much better than a plain round-robin.
    // Balanced routing keeps the natural order and the round-robin.
    int cmax = 0;
    for (int f = 0; f < E; ++f) cmax = max(cmax, s_off[f + 1] - s_off[f]);
    skewed = static_cast<int64_t>(cmax) * E > 2 * static_cast<int64_t>(s_off[E] - s_off[0]);
    for (int e = threadIdx.x; e < E; e += NT) {
      const int c = s_off[e + 1] - s_off[e];
      int r = 0;
      for (int f = 0; f < E; ++f) {
        const int cf = s_off[f + 1] - s_off[f];
        r += (cf > c || (cf == c && f < e)) ? 1 : 0;
      }
      s_tp[skewed ? r : e] = e;
    }
  } else if (warp == 2) {  // tile prefix over experts: ceil(rows / 256)
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int c = e < E ? (s_off[e + 1] - s_off[e] + 2 * BM - 1) / (2 * BM) : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (e < E) s_tp[e] = carry + incl - c;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_tp[E] = carry;
  }
  if (!Tr::kRaggedK && warp == 3) {  // padded offsets: ceil(rows / 128) * 128 per expert
    int carry = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      const int c = e < E ? (s_off[e + 1] - s_off[e] + 127) / 128 * 128 : 0;
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (e < E) s_pad[e] = carry + incl - c;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) s_pad[E] = carry;
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers initialised before any remote arrival
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  const int total = Tr::kRaggedK ? E * p.m_tiles * p.n_tiles : s_tp[E] * p.n_tiles;
  // the it-th tile of this CTA pair (>= total: none left)
  auto tile_at = [&](int it) {
    const int c = (skewed && (it & 1)) ? nclusters - 1 - cluster : cluster;
    return it * nclusters + c;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    // Lane 0 runs the loop alone: no warp collective per stage.
    if (lane == 0) {
      const uint32_t full_cl0 = peer_smem_addr(&full[0], 0);  // CTA 0's full[] (direct mode)
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, arm_par = 0;  // per stage: armed at least once, parity of last arm
      bool ok = true;
      for (int it = 0, tile = tile_at(0); tile < total && ok; tile = tile_at(++it)) {
        const Tile t = decode_tile<MODE>(tile, p, s_tp, s_off, s_pad);
        if constexpr (Tr::kRaggedK) {  // this expert's maps were written by the preceding
          // launch; the thread that issues the copies acquires every map it will use
          if (t.nkb > 0)
            for (int j = 0; j < kMapsPerExpert; ++j) tmap_acquire(p.expert_maps + t.e * kMapsPerExpert + j);
        }
        const int nstage = (t.nkb + HALVES - 1) / HALVES;
        for (int ks = 0; ks < nstage; ++ks) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t *sa = stages + stage * kStageBytes;
          if (rank == 0) {  // both CTAs' bytes
            uint32_t bytes = 2 * kStageBytes;
            if constexpr (!Tr::kRaggedK)
              bytes -= HALVES * (8 - a_boxes(t, 0) - a_boxes(t, 1)) * (32 * BK * 2);
            mbar_arrive_expect_tx(&full[stage], bytes);
          }
          const StageLoad ld{full_cl0 + 8u * stage};
          // a K block past the end (odd count of 64-blocks) loads zero fill or rows
          // that no MMA reads, so every stage carries the same bytes
#pragma unroll
          for (int h = 0; h < HALVES; ++h)
            produce_stage<MODE>(t, ks * HALVES + h, rank, sa + h * kABox, sa + kABytes + h * kBBox, ld,
                                p, &tmA0, &tmA1, &tmB0, &tmB1, &tmA0s, &tmA1s);
          armed |= 1u << stage;
          arm_par = (arm_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      griddep_launch_dependents();  // all loads issued: the next kernel may be launched
      if (*abort_flag && rank == 0) {  // let the pair's copies land before exit
        for (int s = 0; s < STAGES; ++s) {
          if (!((armed >> s) & 1u)) continue;
          for (int i = 0; i < (1 << 22) && !mbar_try_wait(&full[s], (arm_par >> s) & 1u); ++i) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1 && rank == 1) {
    // CTA 1's warp 1 holds the pair's TMEM allocation with CTA 0's warp 1
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (CTA 0)
    // Lane 0 runs the loop alone: no warp collective per stage.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int tile = tile_at(0); tile < total && ok; tile = tile_at(++it)) {
        const Tile t = decode_tile<MODE>(tile, p, s_tp, s_off, s_pad);
        const int buf = it & 1;
        const uint32_t use = (it >> 1) & 1;
        if (!mbar_wait(&tempty[buf], use ^ 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        if (t.nkb == 0) {  // empty expert: both epilogues write zeros
          mbar_arrive(&tfull[buf]);
          mbar_arrive_cluster(peer_smem_addr(&tfull[buf], 1));
          continue;
        }
        const int nstage = (t.nkb + HALVES - 1) / HALVES;
        for (int ks = 0; ks < nstage; ++ks) {
          if (!mbar_wait(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_addr(stages + stage * kStageBytes);
          const uint32_t b_base = a_base + kABytes;
          const int nk16 = (BK / 16) * min(HALVES, t.nkb - ks * HALVES);  // K steps inside K
#pragma unroll
          for (int k16 = 0; k16 < HALVES * (BK / 16); ++k16) {
            if (k16 < nk16) {
              const int h = k16 / (BK / 16), j = k16 % (BK / 16);
              const uint32_t ab = a_base + h * kABox, bb = b_base + h * kBBox;
              const uint64_t adesc = Tr::kAMN ? smem_desc_sw128(ab + j * 2048, kBox, 1024)
                                              : smem_desc_sw128(ab + j * 32, 16, 1024);
              const uint64_t bdesc = Tr::kBMN ? smem_desc_sw128(bb + j * 2048, kBox, 1024)
                                              : smem_desc_sw128(bb + j * 32, 16, 1024);
              tc_mma_f16_pair(d_tmem, adesc, bdesc, Tr::kIdesc, (ks | k16) != 0 ? 1u : 0u);
            }
          }
          tc_commit_pair(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit_pair(&tfull[buf]);
      }
      if (*abort_flag) {  // wait for the pair's MMAs before TMEM is freed
        tc_commit_pair(drain);
        for (int i = 0; i < (1 << 22) && !mbar_try_wait(drain, 0); ++i) {
        }
      }
    }
    __syncwarp();
  } else if (warp < 2 + EW) {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    // column range: warps 2..5 the first, 6..9 the second (a constant 0 with 4 warps)
    const int part = EW == 8 ? (warp - 2) >> 2 : 0;
    const int rit = BM * rank + q * 32 + lane;  // row within the pair's 256-row tile
    const uint32_t tempty0 = peer_smem_addr(&tempty[0], 0);
    const uint32_t tempty1 = peer_smem_addr(&tempty[1], 0);
    // weight quantisation (WQ): the bf16 weight and its codes, [E * wq_rows, wq_ld]
    const int wq_rows = MODE == kFwdGateUp ? p.H : p.I;  // K of the forward GEMM
    const int wq_ld = MODE == kFwdGateUp ? p.I : p.H;
    const SfLayout wq_L{wq_rows, kMxBN};
    const uint16_t *wq_src = p.wsrc[MODE == kFwdGateUp ? rank : 0];
    uint8_t *wq_codes = p.wq[MODE == kFwdGateUp ? rank : 0];
    uint8_t *wq_sf = p.wq_sf[MODE == kFwdGateUp ? rank : 0];
    // The weights for an MXFP8 backward (WQ): of tile i's K blocks (64 weight rows
    // each), the ones of stage ks (128 of K) with ks % (the expert's row tiles)
    // equal to the tile's index among them, so every weight element is quantised
    // once, spread over the expert's tiles.  The epilogue warps share them
    // round-robin in 32-row units and do tile i's after the epilogue of tile
    // i - 1, while tile i's TMA copies bring the same rows into L2, so the
    // weight is read from memory about once.
    auto quant_tile = [&](int i) {
      const int tile = tile_at(i);
      if (tile >= total) return;
      const Tile t = decode_tile<MODE>(tile, p, s_tp, s_off, s_pad);
      const int col0 = MODE == kFwdGateUp ? t.n0 : t.n0 + (BN / 2) * rank;
      if (col0 >= wq_ld) return;
      const int nmt = s_tp[t.e + 1] - s_tp[t.e], mtl = (t.m0 - s_off[t.e]) / (2 * BM);
      int u = 0;
      for (int ks = mtl; ks * HALVES < t.nkb; ks += nmt)
        for (int kb = ks * HALVES; kb < (ks + 1) * HALVES && kb < t.nkb; ++kb)
          for (int q = 0; q < 2; ++q, ++u)
            if ((u + i) % EW == warp - 2)
              quant_weight_rows<MODE == kFwdGateUp ? 4 : 8>(wq_src, t.e * wq_rows + kb * BK + 32 * q, col0,
                                                            wq_ld, wq_codes, wq_sf, wq_L, lane);
    };
    constexpr int kAhead = 1;
    if constexpr (WQ)
      for (int i = 0; i < kAhead; ++i) quant_tile(i);
    int it = 0, gbase = 0;
    for (int tile = tile_at(0); tile < total; tile = tile_at(++it)) {
      const Tile t = decode_tile<MODE>(tile, p, s_tp, s_off, s_pad);
      const int buf = it & 1;
      const uint32_t use = (it >> 1) & 1;
      if (!wait_lane0(&tfull[buf], use, abort_flag)) break;
      __syncwarp();  // every lane reads the accumulator after lane 0 saw it complete
      tc_fence_after();
      const uint32_t tb = tmem_base + buf * BN + (static_cast<uint32_t>(q * 32) << 16);
      uint8_t *stile = epi_tiles + (warp - 2) * kEpiTileBytes;
      if constexpr (MODE == kBwdDA) {
        if (!epilogue_da_ring<Params, BN / 32>(t, tb, rit, q * 32 + lane, p, part, stile, gu_ring,
                                               gu_full, gu_empty, gbase, abort_flag))
          break;
      } else {
        epilogue_tile<MODE>(t, tb, rit, p, part, EW / 4, stile);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(buf ? tempty1 : tempty0);
      if constexpr (WQ) quant_tile(it + kAhead);  // a coming tile's, while its operands stream in
    }
  } else {
    // ------------------------------------------------------------ dA: G/U loader (both CTAs)
    // Walks the tiles in the epilogue's order and loads each tile's G and U,
    // this CTA's 128 rows, in 32-column chunks into the ring (lane 0 alone).
    if (lane == 0) {
      int g = 0;
      uint32_t armed = 0, arm_par = 0;
      bool ok = true;
      for (int it = 0, tile = tile_at(0); tile < total && ok; tile = tile_at(++it)) {
        const Tile t = decode_tile<MODE>(tile, p, s_tp, s_off, s_pad);
        const int nch = min(BN / 32, (p.I - t.n0) / 32);
        for (int c = 0; c < nch; ++c, ++g) {
          const int slot = g % kGuSlots;
          const uint32_t ph = static_cast<uint32_t>(g / kGuSlots) & 1u;
          if (!mbar_wait(&gu_empty[slot], ph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t *dst = gu_ring + slot * kGuChunkBytes;
          mbar_arrive_expect_tx(&gu_full[slot], kGuChunkBytes);
          tma_load_2d(dst, &tmA1, &gu_full[slot], t.n0 + 32 * c, t.m0 + BM * rank);  // G
          tma_load_2d(dst + kGuHalfBytes, &tmB1, &gu_full[slot], t.n0 + 32 * c, t.m0 + BM * rank);  // U
          armed |= 1u << slot;
          arm_par = (arm_par & ~(1u << slot)) | (ph << slot);
        }
      }
      if (*abort_flag) {  // let the copies in flight land before exit
        for (int sl = 0; sl < kGuSlots; ++sl) {
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
  cluster_sync();  // the pair is done with each other's barriers and TMEM
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// Ragged K: per-expert copies of the operand tensor maps whose row extent ends
// at the expert's last row (offsets[e+1]); TMA then zero-fills the rows past it.
struct MapTemplates {
  CUtensorMap m[kMapsPerExpert];
};

__global__ void __launch_bounds__(256) expert_maps_kernel(const __grid_constant__ MapTemplates tm,
                                                          const int32_t *__restrict__ offsets, int E,
                                                          CUtensorMap *out) {
  griddep_wait();  // the previous kernel in the stream has completed
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= E) return;
  const int end = __ldg(offsets + e + 1);
  const uint32_t rows = end > 0 ? static_cast<uint32_t>(end) : 1u;  // an unused map still needs rows >= 1
  for (int j = 0; j < kMapsPerExpert; ++j) {
    const uint4 *src = reinterpret_cast<const uint4 *>(&tm.m[j]);
    CUtensorMap *dst = out + e * kMapsPerExpert + j;
    uint4 *d = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int q = 0; q < 8; ++q) d[q] = src[q];
    tmap_set_global_dim(dst, 1, rows);
  }
  tmap_release();
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// 2-D bf16 tensor map over a row-major [rows, inner] matrix, box {64, box_rows},
// 128-byte swizzle, zero fill out of bounds.
bool make_map(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto fn = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 map over G or U [rows, I]: box {32, 128} (64-byte rows), 64-byte
// swizzle, zero fill out of bounds.
bool make_map_gu(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t rows) {
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

template <int MODE, bool WQ>
cudaError_t launch_kernel(const CUtensorMap &mA0, const CUtensorMap &mA1, const CUtensorMap &mB0,
                          const CUtensorMap &mB1, const CUtensorMap &mA0s, const CUtensorMap &mA1s,
                          const Params &p, int num_sms, cudaStream_t s);

template <int MODE>
cudaError_t launch_mode(const GemmArgs &a, cudaStream_t s) {
  CUtensorMap mA0, mA1, mB0, mB1, mA0s, mA1s;
  Params p{};
  p.M_rows = a.M_rows;
  p.H = a.H;
  p.I = a.I;
  p.E = a.E;
  p.offsets = a.offsets;
  p.o0 = a.o0;
  p.o1 = a.o1;
  p.o2 = a.o2;
  p.o3 = a.o3;
  p.w_row = a.w_row;
  p.aw_t = a.aw_t;
  p.aw_t_sf = a.aw_t_sf;
  p.Mpad = a.Mpad;
  p.g_part = a.g_part;
  p.g_np = 2 * ((a.I + 255) / 256);
  p.status = a.status;
  const uint64_t M = static_cast<uint64_t>(a.M_rows), H = a.H, I = a.I, E = a.E;
  // router modes: a.E is the router's output width, the GEMM sees one expert
  const uint64_t E_out = a.E;
  const bool router = MODE == kRouterFwd || MODE == kRouterDX || MODE == kRouterDW;
  p.E = router ? (MODE == kRouterDW ? (a.r_segments > 0 ? a.r_segments : 1) : 1) : a.E;
  p.of = a.r_out;
  p.n_out = a.E;
  bool ok = true;
  switch (MODE) {
    case kFwdGateUp:
      ok = make_map(&mA0, a.x_perm, H, M, 128) && make_map(&mB0, a.W_gate, I, E * H, 64) &&
           make_map(&mB1, a.W_up, I, E * H, 64) && make_map(&mA0s, a.x_perm, H, M, 32);
      mA1 = mA0;
      mA1s = mA0s;
      p.kdim = a.H;
      p.n_tiles = (a.I + 127) / 128;
      break;
    case kFwdDown:
      ok = make_map(&mA0, a.act, I, M, 128) && make_map(&mB0, a.W_down, H, E * I, 64) &&
           make_map(&mA0s, a.act, I, M, 32);
      mA1 = mA0;
      mA1s = mA0s;
      mB1 = mB0;
      p.kdim = a.I;
      p.n_tiles = (a.H + 255) / 256;
      break;
    case kBwdDA:  // A1, B1: G and U for the epilogue's ring (32 columns x 128 rows)
      ok = make_map(&mA0, a.dy_perm, H, M, 128) && make_map(&mB0, a.W_down, H, E * I, 128) &&
           make_map_gu(&mA1, a.G, I, M) && make_map_gu(&mB1, a.U, I, M) && make_map(&mA0s, a.dy_perm, H, M, 32);
      mA1s = mA0s;
      p.G = a.G;
      p.U = a.U;
      p.kdim = a.H;
      p.n_tiles = (a.I + 255) / 256;
      break;
    case kBwdDX:
      ok = make_map(&mA0, a.dG, I, M, 128) && make_map(&mA1, a.dU, I, M, 128) &&
           make_map(&mB0, a.W_gate, I, E * H, 128) && make_map(&mB1, a.W_up, I, E * H, 128) &&
           make_map(&mA0s, a.dG, I, M, 32) && make_map(&mA1s, a.dU, I, M, 32);
      p.kdim = 2 * a.I;
      p.n_tiles = (a.H + 255) / 256;
      break;
    case kBwdDWDown:
      ok = make_map(&mA0, a.act_w, I, M, 64) && make_map(&mB0, a.dy_perm, H, M, 64);
      mA1 = mA0;
      mB1 = mB0;
      p.m_tiles = (a.I + 2 * BM - 1) / (2 * BM);
      p.n_tiles = (a.H + 255) / 256;
      break;
    case kRouterFwd:  // x [T,H] . W_r [H,E]: one expert, K = H, N = E
      ok = make_map(&mA0, a.r_x, H, M, 128) && make_map(&mB0, a.r_w, E_out, H, 64) &&
           make_map(&mA0s, a.r_x, H, M, 32);
      mA1 = mA0;
      mA1s = mA0s;
      mB1 = mB0;
      p.kdim = a.H;
      p.n_tiles = (a.E + 255) / 256;
      break;
    case kRouterDX:  // bf16(d_logits) [T,E] . W_r^T: K = E (zero-filled to 64s), N = H
      ok = make_map(&mA0, a.r_dlog, E_out, M, 128) && make_map(&mB0, a.r_w, E_out, H, 128) &&
           make_map(&mA0s, a.r_dlog, E_out, M, 32);
      mA1 = mA0;
      mA1s = mA0s;
      mB1 = mB0;
      p.kdim = (a.E + BK - 1) / BK * BK;
      p.n_tiles = (a.H + 255) / 256;
      break;
    case kRouterDW:  // x^T [H,T] . bf16(d_logits) [T,E]: K = T, M = H, N = E
      ok = make_map(&mA0, a.r_x, H, M, 64) && make_map(&mB0, a.r_dlog, E_out, M, 64);
      mA1 = mA0;
      mB1 = mB0;
      p.m_tiles = (a.H + 2 * BM - 1) / (2 * BM);
      p.n_tiles = (a.E + 255) / 256;
      break;
    default:  // kBwdDWGateUp
      ok = make_map(&mA0, a.x_perm, H, M, 64) && make_map(&mB0, a.dG, I, M, 64) &&
           make_map(&mB1, a.dU, I, M, 64);
      mA1 = mA0;
      p.m_tiles = (a.H + 2 * BM - 1) / (2 * BM);
      p.n_tiles = (a.I + 127) / 128;
      break;
  }
  if (!ok) return cudaErrorInvalidValue;
  if constexpr (Traits<MODE>::kRaggedK) {  // whole K blocks: no partial A boxes
    mA0s = mA0;
    mA1s = mA1;
  }
  if constexpr (Traits<MODE>::kRaggedK) {
    if (!a.map_scratch) return cudaErrorInvalidValue;
    MapTemplates tm;
    tm.m[0] = mA0;
    tm.m[1] = mB0;
    tm.m[2] = mB1;
    CUtensorMap *maps = static_cast<CUtensorMap *>(a.map_scratch);
    const cudaError_t e = launch_pdl(expert_maps_kernel, dim3((p.E + 255) / 256), dim3(256), 0, s, 1, tm,
                                     a.offsets, p.E, maps);
    if (e != cudaSuccess) return e;
    p.expert_maps = maps;
  }
  if constexpr (MODE == kFwdGateUp || MODE == kFwdDown) {
    p.wsrc[0] = MODE == kFwdGateUp ? a.W_gate : a.W_down;
    p.wsrc[1] = MODE == kFwdGateUp ? a.W_up : nullptr;
    p.wq[0] = a.wq[0];
    p.wq[1] = a.wq[1];
    p.wq_sf[0] = a.wq_sf[0];
    p.wq_sf[1] = a.wq_sf[1];
    if (a.wq[0]) {  // the variant with weight quantisers
      if (!a.wq_sf[0] || (MODE == kFwdGateUp && (!a.wq[1] || !a.wq_sf[1]))) return cudaErrorInvalidValue;
      return launch_kernel<MODE, true>(mA0, mA1, mB0, mB1, mA0s, mA1s, p, a.num_sms, s);
    }
  }
  return launch_kernel<MODE, false>(mA0, mA1, mB0, mB1, mA0s, mA1s, p, a.num_sms, s);
}

// One launch of a grouped GEMM kernel: clusters of two CTAs, as many pairs as
// fit at once (at most one per two SMs).
template <int MODE, bool WQ>
cudaError_t launch_kernel(const CUtensorMap &mA0, const CUtensorMap &mA1, const CUtensorMap &mB0,
                          const CUtensorMap &mB1, const CUtensorMap &mA0s, const CUtensorMap &mA1s,
                          const Params &p, int num_sms, cudaStream_t s) {
  // once per device: the shared-memory opt-in, and how many CTA pairs fit at once
  static DeviceOnce once;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see launch_pdl
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(threads_of(MODE, WQ));
  cfg.dynamicSmemBytes = smem_bytes(MODE, WQ);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int pair_grid = 0;
  cudaError_t e = once.get(
      [&](int *grid) {
        cudaError_t r = cudaFuncSetAttribute(grouped_gemm_kernel<MODE, WQ>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes(MODE, WQ));
        if (r != cudaSuccess) return r;
        cudaLaunchConfig_t q = cfg;
        q.gridDim = dim3(num_sms & ~1);
        int clusters = 0;
        r = cudaOccupancyMaxActiveClusters(&clusters, grouped_gemm_kernel<MODE, WQ>, &q);
        if (r != cudaSuccess) return r;
        if (clusters < 1) return cudaErrorInvalidConfiguration;
        *grid = 2 * (clusters < num_sms / 2 ? clusters : num_sms / 2);
        return cudaSuccess;
      },
      &pair_grid);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(pair_grid);
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, grouped_gemm_kernel<MODE, WQ>, mA0, mA1, mB0, mB1, mA0s, mA1s, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_grouped_gemm(GemmMode mode, const GemmArgs &a, cudaStream_t s) {
  switch (mode) {
    case kFwdGateUp: return launch_mode<kFwdGateUp>(a, s);
    case kFwdDown: return launch_mode<kFwdDown>(a, s);
    case kBwdDA: return launch_mode<kBwdDA>(a, s);
    case kBwdDX: return launch_mode<kBwdDX>(a, s);
    case kBwdDWDown: return launch_mode<kBwdDWDown>(a, s);
    case kBwdDWGateUp: return launch_mode<kBwdDWGateUp>(a, s);
    case kRouterFwd: return launch_mode<kRouterFwd>(a, s);
    case kRouterDX: return launch_mode<kRouterDX>(a, s);
    case kRouterDW: return launch_mode<kRouterDW>(a, s);
  }
  return cudaErrorInvalidValue;
}

int router_dw_segments(int T, int H, int E) {
  constexpr int kPairs = 76;  // CTA pairs of a 152-SM part
  const int tiles = ((H + 2 * BM - 1) / (2 * BM)) * ((E + 255) / 256);
  int S = kPairs / (tiles > 0 ? tiles : 1);
  S = S < T / 1024 ? S : T / 1024;
  S = S < 32 ? S : 32;
  return S > 1 ? S : 1;
}

const char *gemm_mode_name(GemmMode mode) {
  switch (mode) {
    case kFwdGateUp: return "gemm_gateup_swiglu";
    case kFwdDown: return "gemm_down";
    case kBwdDA: return "gemm_dA_dswiglu";
    case kBwdDX: return "gemm_dX";
    case kBwdDWDown: return "gemm_dW_down";
    case kBwdDWGateUp: return "gemm_dW_gateup";
    case kRouterFwd: return "router_gemm_logits";
    case kRouterDX: return "router_gemm_dx";
    case kRouterDW: return "router_gemm_dW";
  }
  return "?";
}

}  // namespace moe
