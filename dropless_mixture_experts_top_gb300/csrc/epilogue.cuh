// epilogue.cuh -- epilogues of the grouped GEMMs: read one warp's 32 TMEM lanes
// of a 128 x 256 fp32 accumulator and write the layer's bf16 outputs (fused
// SwiGLU for the forward gate/up GEMM, fused dSwiGLU for dA through the G/U
// ring, plain stores for the others, the router projection's fp32 modes).
// epilogue_tile serves both GEMM engines (gemm.cu, and gemm_mx.cu for dX, down
// and the weight gradients; the MXFP8 dA and gate/up epilogues, which also
// quantise, live in gemm_mx.cu).  `P` is any parameter struct with the fields
// used below.
//
// A warp owns 32 rows (one per lane, as tcgen05.ld 32x32b delivers them) and
// walks its columns in 32-column chunks.  Row-major global memory is touched
// through a per-warp 2 KiB shared-memory tile: a lane writes its row's 64
// bytes there, then each instruction moves 8 rows x 64 contiguous bytes
// between the tile and global memory (4 lanes per row), instead of 32 rows x
// 16 bytes.  The tile's 16-byte chunks are XOR-swizzled by row so that both
// access patterns are free of bank conflicts.
#pragma once

#include "common.cuh"
#include "mxfp8.cuh"

namespace moe {

constexpr int kEpiTileBytes = 32 * 32 * 2;  // one warp's 32 x 32 bf16 staging tile

struct Tile {
  int e;        // expert
  int m0;       // first output row of the pair (ragged M: permuted row; ragged K: dW row)
  int row_end;  // ragged M: end of the expert's rows
  int n0;       // first output column
  int nkb;      // K blocks
  int krow0;    // ragged K: expert's first row; ragged M: padded row of m0 (128-aligned segments)
  int kcount;   // ragged K: expert's rows; ragged M: end of the expert's padded segment
};

// Byte offset of row r's 16-byte chunk q (of 4) in a staging tile.
__device__ __forceinline__ uint32_t epi_swz(int r, int q) {
  return static_cast<uint32_t>(r * 64 + ((q ^ ((r >> 1) & 3)) << 4));
}

// The warp's 32 rows x 32 columns, lane = row, to global rows [0, nvalid) at
// g0 (row 0, first column), row stride ld elements.
__device__ __forceinline__ void store_rows32(uint8_t *tile, uint16_t *g0, size_t ld, int nvalid,
                                             const float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
    w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
    w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
    w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
    *reinterpret_cast<uint4 *>(tile + epi_swz(lane, q)) = w;
  }
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 8 * i + (lane >> 2), q = lane & 3;
    const uint4 w = *reinterpret_cast<const uint4 *>(tile + epi_swz(r, q));
    if (r < nvalid) *reinterpret_cast<uint4 *>(g0 + static_cast<size_t>(r) * ld + q * 8) = w;
  }
  __syncwarp();
}

// Coalesced loads of the warp's 32 rows x 32 bf16 columns (rows past nvalid
// read as zero) into registers: issued early, consumed by rows32_to_lanes.
__device__ __forceinline__ void load_rows32(const uint16_t *g0, size_t ld, int nvalid, uint4 (&w)[4]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 8 * i + (lane >> 2), q = lane & 3;
    w[i] = r < nvalid ? __ldg(reinterpret_cast<const uint4 *>(g0 + static_cast<size_t>(r) * ld) + q)
                      : make_uint4(0, 0, 0, 0);
  }
}

// Redistribute loaded rows through the staging tile: lane r gets row r's 32 values.
__device__ __forceinline__ void rows32_to_lanes(uint8_t *tile, const uint4 (&w)[4], float (&v)[32]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = 8 * i + (lane >> 2), q = lane & 3;
    *reinterpret_cast<uint4 *>(tile + epi_swz(r, q)) = w[i];
  }
  __syncwarp();
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 x = *reinterpret_cast<const uint4 *>(tile + epi_swz(lane, q));
    const uint32_t xw[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      v[8 * q + 2 * h] = bf16_lo(xw[h]);
      v[8 * q + 2 * h + 1] = bf16_hi(xw[h]);
    }
  }
  __syncwarp();
}

// The value a bf16 tensor would hold (nearest even), as fp32.
__device__ __forceinline__ float round_bf16(float v) {
  return __uint_as_float(static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v))) << 16);
}

// A warp's 32 x 32 values (lane = row, bf16-exact) quantised down the rows:
// written to the staging tile as bf16, then lane j takes column j's 32 values
// (one 32-token block) and writes its 32 codes at codes + (col0 + j) * ld +
// tok0 and their scale code at sf_byte (its own column's byte).
__device__ __forceinline__ void quant_down_rows32(uint8_t *tile, const float (&v)[32], uint8_t *codes,
                                                  size_t ld, int col0, int tok0, uint8_t *sf_byte) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 w;
    w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
    w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
    w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
    w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
    *reinterpret_cast<uint4 *>(tile + epi_swz(lane, q)) = w;
  }
  __syncwarp();
  float c[32];
  const int qc = lane >> 3, within = (lane & 7) * 2;
#pragma unroll
  for (int i = 0; i < 32; ++i)
    c[i] = __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(
                               tile + epi_swz(i, qc) + within))
                           << 16);
  __syncwarp();  // the tile is rewritten by the next call
  *sf_byte = quant32(c, reinterpret_cast<uint4 *>(codes + static_cast<size_t>(col0 + lane) * ld + tok0));
}

// sigmoid with the approximate (branch-free) reciprocal: within a few fp32 ulp
// of 1 / (1 + e^-z), far below the bf16 rounding of every output it feeds; the
// IEEE division's special-case branch stalled the epilogue warps.
__device__ __forceinline__ float sigmoidf_(float z) { return __fdividef(1.f, 1.f + __expf(-z)); }

__device__ __forceinline__ int clamp_rows(int n) { return n < 0 ? 0 : (n > 32 ? 32 : n); }

// Epilogue of one tile for one warp: 32 rows, and the part-th of nparts column
// ranges (nparts warps share each TMEM lane quarter).  tb: TMEM address of
// this warp's lanes at the accumulator's first column; rit: this lane's row
// within the tile; tile: the warp's staging tile.  NCH: 32-column chunks in
// the tile's unpaired accumulator (8 for 256 columns, 6 for 192); the paired
// modes (gate|up halves) have 4 chunks, each covering both halves.
template <int MODE, class P, int NCH = 8>
__device__ __forceinline__ void epilogue_tile(const Tile &t, uint32_t tb, int rit, const P &p,
                                              int part, int nparts, uint8_t *tile) {
  constexpr int kPairChunks = 4;
  const int cb4 = part * kPairChunks / nparts, ce4 = (part + 1) * kPairChunks / nparts;
  const int cb = part * NCH / nparts, ce = (part + 1) * NCH / nparts;
  const int lane = threadIdx.x & 31;
  uint32_t r0[32], r1[32];
  float v0[32], v1[32], v2[32];
  if constexpr (MODE == kFwdGateUp) {
    const int row = t.m0 + rit, row0 = row - lane;
    const int nvalid = clamp_rows(t.row_end - row0);
    const float w = row < t.row_end ? __ldg(p.w_row + row) : 0.f;
    // for an MXFP8 backward: w * A quantised along tokens -- the warp's 32 rows
    // are one 32-token block of the padded token axis when they start inside
    // the expert's padded segment (rows past its count are zeros)
    const int prow0 = t.krow0 + (rit - lane);
    const bool qtok = p.aw_t != nullptr && prow0 < t.kcount;
    for (int c = cb4; c < ce4; ++c) {
      const int col = t.n0 + 32 * c;
      if (col >= p.I) break;
      tmem_ld32(tb + 32 * c, r0);
      tmem_ld32(tb + 128 + 32 * c, r1);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; i += 2) {  // two columns at a time
        const float g0 = __uint_as_float(r0[i]), g1 = __uint_as_float(r0[i + 1]);
        const float u0 = __uint_as_float(r1[i]), u1 = __uint_as_float(r1[i + 1]);
        const float2 a = f2_get(f2_mul(f2_mul(f2(g0, g1), f2(sigmoidf_(g0), sigmoidf_(g1))), f2(u0, u1)));
        v0[i] = a.x;  // SwiGLU
        v0[i + 1] = a.y;
        v1[i] = g0;
        v1[i + 1] = g1;
        v2[i] = u0;
        v2[i + 1] = u1;
      }
      const size_t off = static_cast<size_t>(row0) * p.I + col;
      store_rows32(tile, p.o0 + off, p.I, nvalid, v0);
      if (p.o1) {  // G, U and w * A are the backward's; a forward that saves nothing skips them
        store_rows32(tile, p.o1 + off, p.I, nvalid, v1);
        store_rows32(tile, p.o2 + off, p.I, nvalid, v2);
      }
      if (p.o3 || qtok) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v0[i] *= w;  // A_w = w * A, the dW_down operand
        if (p.o3) store_rows32(tile, p.o3 + off, p.I, nvalid, v0);
        if (qtok) {  // from the bf16 value the tensor would hold; lane j takes column col + j
          // rows past the count are +0 (0 * A may be -0, whose E4M3 code is not 0)
          const bool valid = row < t.row_end;
#pragma unroll
          for (int i = 0; i < 32; ++i) v1[i] = valid ? round_bf16(v0[i]) : 0.f;
          const int ccol = col + lane;
          const size_t sfb = atom_row_sg<128>(0, ccol, p.Mpad, p.I) + atom_kblock(prow0 >> 5);  // ccol < I: one segment
          quant_down_rows32(tile, v1, p.aw_t, static_cast<size_t>(p.Mpad), col, prow0, p.aw_t_sf + sfb);
        }
      }
    }
  } else if constexpr (MODE == kFwdDown || MODE == kBwdDX) {
    const int row0 = t.m0 + rit - lane;
    const int nvalid = clamp_rows(t.row_end - row0);
    for (int c = cb; c < ce; ++c) {
      const int col = t.n0 + 32 * c;
      if (col >= p.H) break;
      tmem_ld32(tb + 32 * c, r0);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) v0[i] = __uint_as_float(r0[i]);
      store_rows32(tile, p.o0 + static_cast<size_t>(row0) * p.H + col, p.H, nvalid, v0);
    }
  } else if constexpr (MODE == kBwdDWDown) {
    const int i_row0 = t.m0 + rit - lane;
    const int nvalid = clamp_rows(p.I - i_row0);
    for (int c = cb; c < ce; ++c) {
      const int col = t.n0 + 32 * c;
      if (col >= p.H) break;
      if (t.nkb > 0) {
        tmem_ld32(tb + 32 * c, r0);
        tmem_ld_wait();
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) v0[i] = t.nkb > 0 ? __uint_as_float(r0[i]) : 0.f;
      store_rows32(tile, p.o0 + (static_cast<size_t>(t.e) * p.I + i_row0) * p.H + col, p.H, nvalid,
                   v0);
    }
  } else if constexpr (MODE == kRouterFwd || MODE == kRouterDW) {
    // fp32 output [rows, n_out]: logits (rows = tokens, bounded by the segment's
    // end) or dW_r (rows = H, no token ends them; an empty reduction writes 0)
    const int row = t.m0 + rit;
    const bool rv = MODE == kRouterFwd ? row < t.row_end : row < p.H;
    for (int c = cb; c < ce; ++c) {
      const int col = t.n0 + 32 * c;
      if (col >= p.n_out) break;
      if (MODE == kRouterFwd || t.nkb > 0) {
        tmem_ld32(tb + 32 * c, r0);
        tmem_ld_wait();
      }
      if (rv) {  // dW_r split over token segments: segment t.e's partial at t.e * H rows
        const size_t orow = MODE == kRouterDW ? static_cast<size_t>(t.e) * p.H + row : static_cast<size_t>(row);
        float *dst = p.of + orow * p.n_out + col;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (col + 4 * q < p.n_out) {  // n_out is a multiple of 8
            const bool z = MODE == kRouterDW && t.nkb == 0;
            *reinterpret_cast<float4 *>(dst + 4 * q) =
                z ? make_float4(0.f, 0.f, 0.f, 0.f)
                  : make_float4(__uint_as_float(r0[4 * q]), __uint_as_float(r0[4 * q + 1]),
                                __uint_as_float(r0[4 * q + 2]), __uint_as_float(r0[4 * q + 3]));
          }
        }
      }
    }
  } else if constexpr (MODE == kRouterDX) {  // dx [rows, H] bf16 += accumulator
    // K = E is short, so the tile's time is this read-modify-write of dx: the
    // next chunk's rows (other columns) are loaded while this one is processed
    const int row0 = t.m0 + rit - lane;
    const int nvalid = clamp_rows(t.row_end - row0);
    uint16_t *grow = p.o0 + static_cast<size_t>(row0) * p.H;
    uint4 wn[4];
    if (cb < ce && t.n0 + 32 * cb < p.H) load_rows32(grow + t.n0 + 32 * cb, p.H, nvalid, wn);
    for (int c = cb; c < ce; ++c) {
      const int col = t.n0 + 32 * c;
      if (col >= p.H) break;
      uint4 w[4] = {wn[0], wn[1], wn[2], wn[3]};
      uint16_t *g0 = grow + col;
      if (c + 1 < ce && col + 32 < p.H) load_rows32(g0 + 32, p.H, nvalid, wn);
      rows32_to_lanes(tile, w, v1);
      tmem_ld32(tb + 32 * c, r0);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 32; ++i) v0[i] = v1[i] + __uint_as_float(r0[i]);
      store_rows32(tile, g0, p.H, nvalid, v0);
    }
  } else {  // kBwdDWGateUp
    const int h_row0 = t.m0 + rit - lane;
    const int nvalid = clamp_rows(p.H - h_row0);
    for (int c = cb4; c < ce4; ++c) {
      const int col = t.n0 + 32 * c;
      if (col >= p.I) break;
      if (t.nkb > 0) {
        tmem_ld32(tb + 32 * c, r0);
        tmem_ld32(tb + 128 + 32 * c, r1);
        tmem_ld_wait();
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        v0[i] = t.nkb > 0 ? __uint_as_float(r0[i]) : 0.f;
        v1[i] = t.nkb > 0 ? __uint_as_float(r1[i]) : 0.f;
      }
      const size_t off = (static_cast<size_t>(t.e) * p.H + h_row0) * p.I + col;
      store_rows32(tile, p.o0 + off, p.I, nvalid, v0);
      store_rows32(tile, p.o1 + off, p.I, nvalid, v1);
    }
  }
}

// dA's G/U ring (both GEMM engines): a loader warp streams each tile's G and U,
// the CTA's 128 rows, in 32-column chunks (64-byte rows, TMA 64-byte swizzle)
// into kGuSlots slots; the two column halves of epilogue warps take alternate
// chunks, so each half owns one slot.
constexpr int kGuSlots = 2;
constexpr int kGuHalfBytes = 128 * 32 * 2;  // 128 rows x 32 bf16 columns of G (or U): 8 KB
constexpr int kGuChunkBytes = 2 * kGuHalfBytes;

// dA's epilogue for one warp over one tile: its 32 rows, the chunks c of its
// column half (c % 2 == part), G and U taken from the ring that the G/U warp
// fills in chunk order (chunk g of the CTA's sequence sits in slot g %
// kGuSlots; 64-byte rows with the TMA's 64-byte swizzle).  gbase: the CTA's
// running chunk count, advanced past this tile.  With p.g_part set it also
// accumulates the router weight's gradient g_r = <dy_t, Y_r> = <dy_t . W_down^T,
// A_r> over the half's columns (A recomputed from the bf16 G and U, the
// accumulator taken before the router weight) and stores it as partial
// (tile column index, half) of row r.  Returns false if a wait gave up.
template <class P, int NCH>
__device__ __forceinline__ bool epilogue_da_ring(const Tile &t, uint32_t tb, int rit, int rloc,
                                                 const P &p, int part, uint8_t *tile,
                                                 const uint8_t *ring, uint64_t *gu_full,
                                                 uint64_t *gu_empty, int &gbase,
                                                 volatile int *abort_flag) {
  const int lane = threadIdx.x & 31;
  const int row = t.m0 + rit, row0 = row - lane;
  const int nvalid = clamp_rows(t.row_end - row0);
  const float w = row < t.row_end ? __ldg(p.w_row + row) : 0.f;  // dA = w * (dy . W_down^T)
  const size_t rowoff = static_cast<size_t>(row0) * p.I;
  const int nch = min(NCH, (p.I - t.n0) / 32);
  uint32_t r0[32];
  float v1[32], v2[32];
  float gp = 0.f;  // this row's partial router-weight gradient
  bool ok = true;
  for (int c = part; c < nch; c += 2) {
    const int g = gbase + c, slot = g % kGuSlots;
    if (!wait_lane0(&gu_full[slot], static_cast<uint32_t>(g / kGuSlots) & 1u, abort_flag)) {
      ok = false;
      break;
    }
    __syncwarp();  // the other lanes read the chunk after lane 0 saw it land
    const uint8_t *gs = ring + slot * kGuChunkBytes, *us = gs + kGuHalfBytes;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 xg = *reinterpret_cast<const uint4 *>(gs + epi_swz(rloc, q));
      const uint4 xu = *reinterpret_cast<const uint4 *>(us + epi_swz(rloc, q));
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
      const F2 acc = f2(__uint_as_float(r0[i]), __uint_as_float(r0[i + 1]));
      const F2 gg = f2(v1[i], v1[i + 1]), u = f2(v2[i], v2[i + 1]);
      const F2 da = f2_mul(w2, acc);
      const F2 sg = f2(sigmoidf_(v1[i]), sigmoidf_(v1[i + 1]));
      const F2 silu = f2_mul(gg, sg);
      const float2 su = f2_get(f2_mul(silu, u));
      gp = fmaf(__uint_as_float(r0[i]), su.x, gp);  // <dy . W_down^T, A>, in column order
      gp = fmaf(__uint_as_float(r0[i + 1]), su.y, gp);
      const float2 dg = f2_get(f2_mul(f2_mul(f2_mul(da, u), sg), f2_fma(gg, f2_sub(one, sg), one)));
      const float2 du = f2_get(f2_mul(da, silu));  // dU = dA * silu(G)
      v2[i] = dg.x;
      v2[i + 1] = dg.y;
      v1[i] = du.x;
      v1[i + 1] = du.y;
    }
    store_rows32(tile, p.o0 + rowoff + col, p.I, nvalid, v2);
    store_rows32(tile, p.o1 + rowoff + col, p.I, nvalid, v1);
  }
  if (ok && p.g_part && row < t.row_end)
    p.g_part[static_cast<size_t>(row) * p.g_np + (t.n0 >> 8) * 2 + part] = gp;
  gbase += nch;
  return ok;
}

}  // namespace moe
